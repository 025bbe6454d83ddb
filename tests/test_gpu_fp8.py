"""fp8 (E4M3) KV cache on the GPU, through the C ABI, against the oracle:
the quantizing append and the block copy bit for bit, attention over E4M3
pools within the attention tolerance. Pool rows no sequence may read hold the
E4M3 NaN code, so a read outside a sequence's tokens fails the comparison."""

import math

import numpy as np
import pytest

import oracle
import synthetic
from tests.gpu_helpers import assert_close_attention, used_rows_mask

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

NAN8 = np.uint8(0x7F)


@pytest.fixture(scope="module")
def pa(libpa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return libpa


def d(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _scales(rng, hkv):
    return (rng.uniform(0.002, 0.02, hkv).astype(np.float32),
            rng.uniform(0.002, 0.02, hkv).astype(np.float32))


def _fp8_case(seed, S, Hq, Hkv, D, BS, lens, nb_extra=3):
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
    kp = synthetic.fp8_codes(rng, (nb, BS, Hkv, D))
    vp = synthetic.fp8_codes(rng, (nb, BS, Hkv, D))
    keep = used_rows_mask(table, lens, nb, BS)
    kp[~keep] = NAN8
    vp[~keep] = NAN8
    ks, vs = _scales(rng, Hkv)
    return q, kp, vp, ks, vs, table


def _attend(pa, q, kp, vp, ks, vs, table, lens, scale, partition=0):
    out = pa.pa_decode_attention_fp8(d(q), d(kp), d(vp), d(ks), d(vs), d(table.astype(np.int32)),
                                     d(np.asarray(lens, np.int32)), scale,
                                     partition_tokens=partition)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_append_fp8_bit_exact(pa):
    rng = np.random.default_rng(21)
    NB, BS, H, D = 9, 16, 4, 128
    kp = synthetic.fp8_codes(rng, (NB, BS, H, D))
    vp = synthetic.fp8_codes(rng, (NB, BS, H, D))
    T = 12
    kn = (rng.standard_normal((T, H, D)) * 3).astype(np.float16)
    vn = (rng.standard_normal((T, H, D)) * 3).astype(np.float16)
    # saturation, subnormal and zero codes must come out exactly too
    kn[0, 0, :8] = np.array([60000, -60000, 1e-4, -1e-4, 0, -0.0, 5e-3, 7.0], np.float16)
    vn[1, 2, :4] = np.array([-30000, 2e-5, 0, 3.5], np.float16)
    ks, vs = _scales(rng, H)
    slots = np.array([0, 17, 35, -1, 143, 100, 5, 63, 64, 80, -1, 15], np.int32)
    dk, dv = d(kp), d(vp)
    pa.pa_append_kv_fp8(d(kn), d(vn), dk, dv, d(slots), d(ks), d(vs))
    torch.cuda.synchronize()
    ek, ev = oracle.append_kv_fp8(kp, vp, kn, vn, slots, ks, vs)
    assert np.array_equal(dk.cpu().numpy(), ek)
    assert np.array_equal(dv.cpu().numpy(), ev)
    assert pa.pa_device_error() == 0


def test_copy_blocks_fp8_bit_exact(pa):
    rng = np.random.default_rng(22)
    NB, BS, H, D = 8, 16, 2, 128
    kp = rng.integers(0, 256, (NB, BS, H, D), dtype=np.uint8)
    vp = rng.integers(0, 256, (NB, BS, H, D), dtype=np.uint8)
    pairs = np.array([[1, 4], [6, 0], [2, 7]], np.int32)
    dk, dv = d(kp), d(vp)
    pa.pa_copy_blocks_fp8(dk, dv, d(pairs))
    torch.cuda.synchronize()
    ek, ev = oracle.copy_blocks(kp, vp, pairs)
    assert np.array_equal(dk.cpu().numpy(), ek)
    assert np.array_equal(dv.cpu().numpy(), ev)


@pytest.mark.parametrize("BS", [16, 32])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_fp8_shape_matrix(pa, BS, G):
    Hkv = 2
    lens = [1, BS - 1, BS, BS + 1, 255, 256, 257, 700]
    q, kp, vp, ks, vs, table = _fp8_case(BS * 10 + G, len(lens), G * Hkv, Hkv, 128, BS, lens)
    scale = np.float32(1 / math.sqrt(128))
    got = _attend(pa, q, kp, vp, ks, vs, table, lens, scale)
    exp = oracle.decode_attention_fp8(q, kp, vp, ks, vs, table, lens, scale)
    assert_close_attention(got, exp, f"fp8 BS{BS} G{G}")
    assert pa.pa_device_error() == 0


@pytest.mark.parametrize("partition", [16, 48, 256])
def test_fp8_partitions(pa, partition):
    lens = [1, 300, 1000, 4097]
    q, kp, vp, ks, vs, table = _fp8_case(31, 4, 16, 4, 128, 16, lens)
    got = _attend(pa, q, kp, vp, ks, vs, table, lens, np.float32(0.088), partition)
    exp = oracle.decode_attention_fp8(q, kp, vp, ks, vs, table, lens, np.float32(0.088))
    assert_close_attention(got, exp, f"fp8 partition {partition}")


def test_fp8_zero_length(pa):
    lens = [0, 5, 0, 40]
    q, kp, vp, ks, vs, table = _fp8_case(32, 4, 8, 2, 128, 16, [1, 5, 1, 40])
    got = _attend(pa, q, kp, vp, ks, vs, table, lens, np.float32(0.1))
    assert not got[0].any() and not got[2].any()
    exp = oracle.decode_attention_fp8(q, kp, vp, ks, vs, table, lens, np.float32(0.1))
    assert_close_attention(got, exp, "fp8 zero length")


@pytest.mark.parametrize("every_code", [False, True])
def test_fp8_gqa_batch_full_size_sampled(pa, every_code):
    """The 64-sequence GQA batch (lengths U[128, 2048], 32q/8kv, D=128,
    BS=16) over an E4M3 cache, in the launch configuration the benchmark
    uses; every head of sampled sequences checked against the oracle. The
    cache's codes are those of a scaled N(0,1) tensor, or every finite code
    equally often (zeros, subnormals, every exponent field, +-448)."""
    b = synthetic.config2_gqa_batch()
    c = synthetic.fp8_cache(b, every_code=every_code)
    ref = oracle.decode_step(b, compute_attention=False)
    keep = used_rows_mask(ref.block_table, ref.seq_lens, b.num_blocks, b.block_size)
    kp, vp = c.k_pool.copy(), c.v_pool.copy()
    kp[~keep] = NAN8
    vp[~keep] = NAN8
    got = _attend(pa, b.q, kp, vp, c.k_scale, c.v_scale, ref.block_table, ref.seq_lens, b.scale)
    seqs = [0, 17, 40, 63]
    exp = oracle.decode_attention_fp8(b.q, kp, vp, c.k_scale, c.v_scale, ref.block_table,
                                      ref.seq_lens, b.scale, seqs=seqs)
    assert_close_attention(got[seqs], exp[seqs], "fp8 gqa batch")
    assert np.isfinite(got).all()


def test_fp8_append_then_attend(pa):
    """One decode step on an E4M3 cache: quantizing append of the new token,
    then attention over every cached token including it."""
    rng = np.random.default_rng(40)
    lens_before = [30, 15, 200]
    S, Hq, Hkv, D, BS = 3, 8, 2, 128, 16
    lens = [L + 1 for L in lens_before]
    q, kp, vp, ks, vs, table = _fp8_case(41, S, Hq, Hkv, D, BS, lens)
    slots = np.array([int(table[i, L // BS]) * BS + L % BS for i, L in enumerate(lens_before)],
                     np.int32)
    kn = rng.standard_normal((S, Hkv, D)).astype(np.float16)
    vn = rng.standard_normal((S, Hkv, D)).astype(np.float16)
    dk, dv = d(kp), d(vp)
    pa.pa_append_kv_fp8(d(kn), d(vn), dk, dv, d(slots), d(ks), d(vs))
    out = pa.pa_decode_attention_fp8(d(q), dk, dv, d(ks), d(vs), d(table), d(np.asarray(lens, np.int32)),
                                     np.float32(0.09))
    torch.cuda.synchronize()
    ek, ev = oracle.append_kv_fp8(kp, vp, kn, vn, slots, ks, vs)
    assert np.array_equal(dk.cpu().numpy(), ek) and np.array_equal(dv.cpu().numpy(), ev)
    exp = oracle.decode_attention_fp8(q, ek, ev, ks, vs, table, lens, np.float32(0.09))
    assert_close_attention(out.cpu().numpy(), exp, "fp8 step")


@pytest.mark.parametrize("D,BS", [(64, 16), (128, 8)])
def test_fp8_unsupported_shapes_are_refused(pa, D, BS):
    from paged_kv_cache_40_gb300 import PaError
    lens = [20]
    q, kp, vp, ks, vs, table = _fp8_case(50, 1, 2, 2, D, BS, lens)
    with pytest.raises(PaError):
        _attend(pa, q, kp, vp, ks, vs, table, lens, np.float32(0.1))


# ---------------------------------------------------- every finite E4M3 code --
def _every_code_case(seed, lens, G, Hkv, BS):
    """Pools whose attended rows hold every finite E4M3 code (each equally
    often, seeded order) and whose other rows hold the NaN code."""
    rng = np.random.default_rng(seed)
    S, D = len(lens), 128
    mb = max(1, max(-(-L // BS) for L in lens))
    nb = sum(-(-L // BS) for L in lens) + 3
    perm = rng.permutation(nb)
    table = -np.ones((S, mb), np.int32)
    pos = 0
    for i, L in enumerate(lens):
        n = -(-L // BS)
        table[i, :n] = perm[pos:pos + n]
        pos += n
    keep = used_rows_mask(table, lens, nb, BS)
    kp = np.full((nb, BS, Hkv, D), NAN8, np.uint8)
    vp = np.full((nb, BS, Hkv, D), NAN8, np.uint8)
    rows = int(keep.sum())
    kp[keep] = synthetic.fp8_codes_every_finite(rng, (rows, Hkv, D))
    vp[keep] = synthetic.fp8_codes_every_finite(rng, (rows, Hkv, D))
    finite = set(synthetic.fp8_finite_codes().tolist())
    assert set(np.unique(kp[keep]).tolist()) == finite
    assert set(np.unique(vp[keep]).tolist()) == finite
    q = rng.standard_normal((S, G * Hkv, D)).astype(np.float16)
    ks, vs = _scales(rng, Hkv)
    return q, kp, vp, ks, vs, table


@pytest.mark.parametrize("layout", ["pools", "records"])
@pytest.mark.parametrize("BS", [16, 32])
@pytest.mark.parametrize("G", [1, 4, 8])
def test_fp8_every_finite_code(pa, layout, BS, G):
    """Attention over E4M3 pools holding every finite code (zero and -0,
    +-subnormals, exponent fields 1..15, the saturation value +-448), in two
    pools and in the one-pool record layout, against the oracle's attention
    of the decoded values."""
    lens = [1, BS - 1, BS, BS + 1, 300, 777]
    Hkv = 2
    q, kp, vp, ks, vs, table = _every_code_case(600 + 10 * BS + G, lens, G, Hkv, BS)
    scale = np.float32(1 / math.sqrt(128))
    if layout == "pools":
        got = _attend(pa, q, kp, vp, ks, vs, table, lens, scale)
        exp = oracle.decode_attention_fp8(q, kp, vp, ks, vs, table, lens, scale)
    else:
        recs = oracle.make_kv_pool(kp, vp)
        raw = recs.view(np.uint8).reshape(len(recs), 2, BS, Hkv, 128)
        kv = d(raw)
        k, v = pa.kv_views(kv)
        out = pa.pa_decode_attention_fp8(d(q), k, v, d(ks), d(vs), d(table),
                                         d(np.asarray(lens, np.int32)), scale)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        exp = oracle.decode_attention_interleaved_fp8(q, recs, ks, vs, table, lens, scale)
    assert np.isfinite(got).all()
    assert_close_attention(got, exp, f"fp8 every code {layout} BS{BS} G{G}")
    assert pa.pa_device_error() == 0
