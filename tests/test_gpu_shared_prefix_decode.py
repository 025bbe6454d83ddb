"""pa_decode_attention_shared_prefix on the GPU (through the C ABI) against the
fp64 oracle's plain attention: sequences that share their first P physical
blocks, with private suffixes of every length class. Rows no sequence may read
are NaN-poisoned."""

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


def d(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _case(seed, S, Hq, Hkv, BS, P, suffix_lens, D=128, extra=4, mb=None):
    """P shared blocks, then per-sequence private blocks for its suffix; the
    table is P + the longest suffix's blocks + 1 wide unless `mb` is given."""
    rng = np.random.default_rng(seed)
    lens = [P * BS + s for s in suffix_lens]
    priv = [-(-s // BS) for s in suffix_lens]
    nb = P + sum(priv) + extra
    perm = rng.permutation(nb).astype(np.int32)
    prefix = perm[:P]
    mb = P + max(priv) + 1 if mb is None else mb
    table = -np.ones((S, mb), np.int32)
    pos = P
    for i in range(S):
        table[i, :P] = prefix
        table[i, P:P + priv[i]] = perm[pos:pos + priv[i]]
        pos += priv[i]
    q = rng.standard_normal((S, Hq, D)).astype(np.float16)
    kp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    vp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    kp, vp = poison_unread_rows(kp, vp, table, lens, BS)
    return q, kp, vp, prefix, table, np.asarray(lens, np.int32)


def _run(pa, q, kp, vp, prefix, table, lens, scale):
    out = pa.pa_decode_attention_shared_prefix(d(q), d(kp), d(vp), d(prefix), d(table), d(lens),
                                               scale)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("BS", [16, 32])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_shared_prefix_matrix(pa, BS, G):
    Hkv = 2
    suffix = [0, 1, BS - 1, BS, 3 * BS + 5, 200, 7]
    q, kp, vp, prefix, table, lens = _case(BS * 10 + G, len(suffix), G * Hkv, Hkv, BS, 5, suffix)
    scale = np.float32(1 / math.sqrt(128))
    got = _run(pa, q, kp, vp, prefix, table, lens, scale)
    exp = oracle.decode_attention(q, kp, vp, table, lens, scale)
    assert_close_attention(got, exp, f"shared prefix BS{BS} G{G}")
    assert pa.pa_device_error() == 0


def test_shared_prefix_many_rows_and_chunks(pa):
    """300 sequences (19 row tiles of 64 (sequence, head) rows per KV head)
    over a 96-block prefix split into chunks."""
    rng = np.random.default_rng(3)
    suffix = rng.integers(0, 80, 300).tolist()
    q, kp, vp, prefix, table, lens = _case(4, 300, 32, 8, 16, 96, suffix)
    got = _run(pa, q, kp, vp, prefix, table, lens, np.float32(0.088))
    seqs = [0, 1, 63, 64, 150, 299]
    exp = oracle.decode_attention(q, kp, vp, table, lens, np.float32(0.088), seqs=seqs)
    assert_close_attention(got[seqs], exp[seqs], "many rows")
    assert np.isfinite(got).all()


def test_shared_prefix_first_step_of_prefix_workload(pa):
    """The shared-prefix workload's first decode step (128 sequences forked
    from one 2040-token prefix, 32q/8kv): tables from the native block
    manager after the copy-on-write step; the 127 full prefix blocks are the
    shared prefix."""
    w = synthetic.config4_shared_prefix()
    a = pa.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    a.add_seq(0, w.prefix_len)
    for c in range(1, w.num_seqs):
        a.fork(0, c)
    active = list(range(w.num_seqs))
    a.append_slots(active)
    mb = -(-(w.prefix_len + 1) // w.block_size)
    table, lens = a.build_tables(active, mb)
    P = w.prefix_len // w.block_size
    prefix = table[0, :P].copy()
    assert (table[:, :P] == prefix).all()
    q = w.step_inputs(0, w.num_seqs)[0]
    got = _run(pa, q, w.k_pool, w.v_pool, prefix, table, lens, w.scale)
    seqs = [0, 5, 64, 127]
    exp = oracle.decode_attention(q, w.k_pool, w.v_pool, table, lens, w.scale, seqs=seqs)
    assert_close_attention(got[seqs], exp[seqs], "prefix workload first step")


def test_zero_prefix_blocks_is_plain_decode(pa):
    q, kp, vp, prefix, table, lens = _case(8, 3, 8, 2, 16, 0, [5, 40, 300])
    got = _run(pa, q, kp, vp, np.zeros(0, np.int32), table, lens, np.float32(0.1))
    exp = oracle.decode_attention(q, kp, vp, table, lens, np.float32(0.1))
    assert_close_attention(got, exp, "P = 0")


def test_sequence_shorter_than_prefix_is_reported(pa):
    q, kp, vp, prefix, table, lens = _case(9, 2, 8, 2, 16, 4, [3, 3])
    lens = lens.copy()
    lens[1] = 20                                   # 4 prefix blocks hold 64 tokens
    _run(pa, q, kp, vp, prefix, table, lens, np.float32(0.1))
    with pytest.raises(pa.PaError) as e:
        pa.pa_device_error()
    assert e.value.flags & pa.PA_DEVERR_BAD_LEN


# ------------------------------------------------ short suffixes: one launch --
# A table at most 32 tokens wider than the prefix means every suffix is that
# short: the call then runs as one launch whose clusters (the prefix chunks of
# a row tile and KV head) merge their partials on chip and attend the
# suffixes themselves. Cluster sizes 8, 4, 2 and 1 come from the prefix
# length and the grid; chunks past a short prefix are empty.
@pytest.mark.parametrize("BS", [16, 32])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("P", [1, 2, 5, 9])
def test_short_suffix_one_launch_matrix(pa, BS, G, P):
    Hkv = 2
    suffix = [0, 1, 7, BS - 1, BS, 32, 31, 2, 0, 17, 32]
    q, kp, vp, prefix, table, lens = _case(1000 + 100 * P + BS + G, len(suffix), G * Hkv, Hkv,
                                           BS, P, suffix, mb=P + 32 // BS)
    scale = np.float32(1 / math.sqrt(128))
    got = _run(pa, q, kp, vp, prefix, table, lens, scale)
    exp = oracle.decode_attention(q, kp, vp, table, lens, scale)
    assert_close_attention(got, exp, f"short suffix BS{BS} G{G} P{P}")
    assert pa.pa_device_error() == 0


@pytest.mark.parametrize("S,G,Hkv", [(128, 4, 8), (300, 4, 8), (40, 8, 8), (3, 1, 1)])
def test_short_suffix_one_launch_grids(pa, S, G, Hkv):
    """Row tiles x KV heads x cluster sizes across the grid's range: the
    prefix workload's shape (4 row tiles, clusters of 4), 10 row tiles (no
    cluster), one row tile of 8 heads, a single row."""
    rng = np.random.default_rng(S)
    suffix = rng.integers(0, 17, S).tolist()
    P = 40
    q, kp, vp, prefix, table, lens = _case(7 + S, S, G * Hkv, Hkv, 16, P, suffix, mb=P + 1)
    got = _run(pa, q, kp, vp, prefix, table, lens, np.float32(0.088))
    seqs = sorted({0, 1, S // 2, S - 1})
    exp = oracle.decode_attention(q, kp, vp, table, lens, np.float32(0.088), seqs=seqs)
    assert_close_attention(got[seqs], exp[seqs], f"short suffix S{S} G{G} Hkv{Hkv}")
    assert np.isfinite(got).all()
    assert pa.pa_device_error() == 0


def test_short_suffix_bad_length_and_block_are_reported(pa):
    q, kp, vp, prefix, table, lens = _case(11, 4, 8, 2, 16, 6, [3, 9, 16, 0], mb=8)
    lens = lens.copy()
    lens[3] = 6 * 16 - 5                           # shorter than the prefix
    _run(pa, q, kp, vp, prefix, table, lens, np.float32(0.1))
    with pytest.raises(pa.PaError) as e:
        pa.pa_device_error()
    assert e.value.flags & pa.PA_DEVERR_BAD_LEN
    table = table.copy()
    table[1, 6] = 10_000_000                       # a suffix block outside the pool
    lens[3] = 6 * 16
    _run(pa, q, kp, vp, prefix, table, lens, np.float32(0.1))
    with pytest.raises(pa.PaError) as e:
        pa.pa_device_error()
    assert e.value.flags & pa.PA_DEVERR_BAD_BLOCK


# ---------------------------------- short suffixes on the tensor cores --
# In the one-launch mode the CTA that finishes a slice of a tile's rows also
# attends the suffixes of that slice's sequences, as extra 128-token
# sub-chunks: W = (table width - P) * BS tokens per sequence, 128 / W
# sequences per sub-chunk, each row masked to its own sequence's tokens; V
# rows past a length are cleared before the P V MMAs (the poisoned rows here
# would otherwise reach the output as 0 * NaN).
@pytest.mark.parametrize("scale", [0.088, -0.07, 0.6])
def test_two_suffix_subchunks_and_an_empty_chunk(pa, scale):
    """64 sequences, G = 2: one row tile in clusters of 4 chunks over a
    5-block prefix (the last chunk holds no prefix block), 16 sequences per
    slice with 16 suffix tokens each = two suffix sub-chunks per CTA; the
    last CTA's rows have only suffix sub-chunks. At scale 0.6 the running
    max often moves by more than 2^8, so O is rescaled in tensor memory."""
    rng = np.random.default_rng(21)
    suffix = rng.integers(0, 17, 64).tolist()
    suffix[:4] = [0, 16, 1, 15]
    suffix[-3:] = [0, 16, 3]
    q, kp, vp, prefix, table, lens = _case(31, 64, 4, 2, 16, 5, suffix, mb=6)
    got = _run(pa, q, kp, vp, prefix, table, lens, np.float32(scale))
    exp = oracle.decode_attention(q, kp, vp, table, lens, np.float32(scale))
    assert_close_attention(got, exp, f"two suffix sub-chunks, scale {scale}")
    assert pa.pa_device_error() == 0


def test_suffix_width_32_in_two_subchunks(pa):
    """128 sequences, 32 q / 8 kv heads, a 40-block prefix and a table two
    blocks wider: 8 sequences per slice x 32 suffix tokens = two sub-chunks."""
    rng = np.random.default_rng(22)
    suffix = rng.integers(0, 33, 128).tolist()
    suffix[:5] = [0, 32, 16, 17, 31]
    q, kp, vp, prefix, table, lens = _case(32, 128, 32, 8, 16, 40, suffix, mb=42)
    got = _run(pa, q, kp, vp, prefix, table, lens, np.float32(0.088))
    seqs = [0, 1, 2, 3, 4, 63, 64, 127]
    exp = oracle.decode_attention(q, kp, vp, table, lens, np.float32(0.088), seqs=seqs)
    assert_close_attention(got[seqs], exp[seqs], "suffix width 32")
    assert np.isfinite(got).all()
    assert pa.pa_device_error() == 0


def test_zero_scale_gives_uniform_weights(pa):
    """scale 0: every token of a sequence weighs the same (the call takes the
    two-kernel path for it)."""
    suffix = [0, 1, 9, 16, 5]
    q, kp, vp, prefix, table, lens = _case(33, 5, 8, 2, 16, 6, suffix, mb=7)
    got = _run(pa, q, kp, vp, prefix, table, lens, np.float32(0.0))
    exp = oracle.decode_attention(q, kp, vp, table, lens, np.float32(0.0))
    assert_close_attention(got, exp, "scale 0")
    assert pa.pa_device_error() == 0
