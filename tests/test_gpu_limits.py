"""Decode attention at the limits of what the library serves, on the GPU
against the oracle: the largest batch (16384 sequences, the prefix sum over
all of them in shared memory), and the degenerate batch in which no sequence
has a token. Unread pool rows are NaN-poisoned."""

import numpy as np
import pytest

import oracle
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


def _batch(seed, lens, Hq, Hkv, D, BS):
    rng = np.random.default_rng(seed)
    S = len(lens)
    mb = max(1, max(-(-int(L) // BS) for L in lens))
    nb = sum(-(-int(L) // BS) for L in lens) + 3
    perm = rng.permutation(nb).astype(np.int32)
    table = -np.ones((S, mb), np.int32)
    pos = 0
    for i, L in enumerate(lens):
        n = -(-int(L) // BS)
        table[i, :n] = perm[pos:pos + n]
        pos += n
    q = rng.standard_normal((S, Hq, D)).astype(np.float16)
    kp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    vp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    kp, vp = poison_unread_rows(kp, vp, table, lens, BS)
    return q, kp, vp, table


def test_largest_batch_16384_sequences(pa):
    rng = np.random.default_rng(77)
    S = 16384
    lens = rng.integers(0, 41, S).astype(np.int32)
    lens[[5, 16383]] = 0
    lens[[0, 8191]] = 40
    q, kp, vp, table = _batch(78, lens, 8, 2, 64, 16)
    out = pa.pa_decode_attention(d(q), d(kp), d(vp), d(table), d(lens), np.float32(0.125))
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert pa.pa_device_error() == 0
    assert np.isfinite(got).all()
    assert not got[5].any() and not got[16383].any()
    seqs = [0, 1, 2, 777, 8191, 8192, 12000, 16382] + rng.integers(0, S, 8).tolist()
    exp = oracle.decode_attention(q, kp, vp, table, lens, np.float32(0.125), seqs=seqs)
    assert_close_attention(got[seqs], exp[seqs], "16384 sequences")


def test_batch_with_no_tokens_at_all(pa):
    q, kp, vp, table = _batch(79, [1, 1, 1, 1, 1], 8, 2, 128, 16)
    lens = np.zeros(5, np.int32)
    out = torch.full(q.shape, 7.0, dtype=torch.float16, device="cuda")
    pa.pa_decode_attention(d(q), d(kp), d(vp), d(table), d(lens), 0.1, out=out)
    torch.cuda.synchronize()
    assert not out.any()
    assert pa.pa_device_error() == 0
